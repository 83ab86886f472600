// qmv_mtile.cu -- M-column tiles on the bulk-copy pipeline (M >= 2 token
// columns, K a multiple of 256).
//
// What they compute ("raw-metal-loop-playbook", prefill-regimes table: keep
// each output scalar's K-dot in the single-token accumulation order and stage
// the weights across the M columns): every column is bit-identical to the
// M = 1 pipeline's result for that column, in the exact form (the oracle's
// order) and in the fast mode's folded-offset form (see qmv_decode.cuh) --
// the same per-block chains, block finish and serial fold over the blocks.
//
// Layout of the work:
//   * a segment's activation table depends on the activations only, not on
//     the weight rows, so a small kernel first builds every (column chunk,
//     512-code segment) table once per call, with its block sums, into the
//     caller's workspace (8960 bytes each for 4 columns, 17408 for 8; a few
//     hundred KB that stay in L2);
//   * a tile is R = 32*U weight rows x MC = 4 or 8 token columns over the
//     whole K (a cost model picks U and MC; with 8 columns each code's mask
//     serves twice the paired FMAs, and two ring stages fit); a persistent
//     CTA (one per SM) walks its tiles, each in segments of 512 codes;
//   * the copy warp brings, per segment, the tile's packed codes (one or more
//     128-byte-swizzled boxes of R rows x 128 bytes), its group-32 scales and
//     the segment's prebuilt table into a ring of stages;
//   * each 64-code item of the segment goes to one compute warp (two for
//     128-row, 4-column tiles, each taking half the rows): lane l holds rows
//     l + 32u,
//     decodes each code once and runs the paired-FMA chains of the MC columns
//     (one 16-byte shared-memory broadcast serves two columns of its rows);
//     the block results go to one of two fold buffers (one 16-byte store per
//     row), so the compute warps only decode and FMA;
//   * the fold warps (four, or two beside sixteen compute warps), one segment
//     behind, add the block results in block order: each thread owns some
//     rows' (row, column) accumulators, and stores them after the tile's last
//     segment.
// With the fused residual-add + RMSNorm prologue, the table kernel forms
// each of its columns' h = fp16(x + r), the sum of squares in the oracle's
// order and inv, then the normalised fp16 activations y = fp16((h*inv)*gamma)
// of its segment, from which it builds the table, and stores that segment of
// h to h_out: once per column and segment instead of once per row tile, and
// y is what the fused definition feeds the matvec.
// The roles meet only on mbarriers (stage full/empty, fold buffer
// full/empty), so a slow warp delays the others by its lag, not by a
// CTA-wide barrier per segment.  Every wait is bounded; a wait that runs out
// records an error code in this file's device error word and the CTA winds
// down.
#include <cuda.h>

#include "qmv_pipe.cuh"
#include "qmv_prologue.cuh"

namespace qmv {

__device__ int g_mt_error = 0;

namespace {

using namespace pipe;

constexpr int MT_NSMAX = 3;                  // ring stages (at most)
constexpr int MT_KS = 512;                   // codes per segment
constexpr int MT_ITEMS = MT_KS / 64;         // 64-code items per segment (one per compute warp)
constexpr int MT_BLOCKS = MT_KS / 32;        // 32-code blocks per segment
constexpr int MT_HDR = 1024;                 // barriers, flags
constexpr int ERR_MT_TIMEOUT = 32;

// One segment's table record for MC token columns, as the table kernel
// writes it to the workspace and the copy warp brings it into a stage: per
// item 4 octets of 8 steps, a step MC fp32 pairs (the columns side by side),
// each octet padded by 16 bytes, then the block sums [block][MC] (fast mode).
template <int MC>
struct MtRec {
  static constexpr int OCT = 8 * MC + 2;                 // u64 per octet
  static constexpr int TITEM = 4 * OCT;                  // u64 per item
  static constexpr int TAB = MT_ITEMS * TITEM * 8;       // table bytes
  static constexpr int YSUM = MT_BLOCKS * MC * 4;        // block-sum bytes
  static constexpr int TBLK = TAB + YSUM;                // 8960 (MC 4) or 17408 (MC 8) bytes
  static_assert(TBLK % 256 == 0, "records start 256-byte aligned in the workspace; bulk copies move 16-byte multiples");
};
constexpr int MT_TB_THREADS = 32;                        // threads of the table kernel per column

// Shared-memory layout of one kernel variant (offsets from a 1024-byte
// aligned base; the copies with 128-byte swizzle need 1024-byte aligned
// boxes).
template <int BITS, int U, int MC_>
struct MtLayout {
  static constexpr int MC = MC_;                           // token columns per tile (4 or 8)
  static constexpr int R = 32 * U;                         // rows per tile
  static constexpr int NS = (MC == 8) ? 2 : 3;             // ring stages (what fits)
  static constexpr int TBLK = MtRec<MC>::TBLK;
  // 128-row tiles of 4 columns split each item's rows over two compute warps
  // (four per scheduler: more warps to hide the paired FMAs' and loads'
  // latencies); other tiles keep one warp per item (their FMA chains are
  // long enough, or their rows are few)
  static constexpr int CWI = (U >= 4 && MC == 4) ? 2 : 1;  // compute warps per item (row halves)
  static constexpr int UW = U / CWI;                       // rows per lane of a compute warp
  static constexpr int CW = MT_ITEMS * CWI;                // compute warps
  static constexpr int TW = (CWI == 2) ? 2 : 4;            // fold warps (within the register file)
  static constexpr int THREADS = 32 * (CW + TW + 1);       // + fold warps + the copy warp
  static constexpr int NBOX = BITS / 2;                    // 128-byte code boxes per row per segment
  static constexpr int BOX = R * 128;
  static constexpr int SC_OFF = NBOX * BOX;                // scales: [R][16] fp16
  static constexpr int TBL_OFF = SC_OFF + R * 32;          // the segment's table record
  static constexpr int STAGE = (TBL_OFF + TBLK + 1023) / 1024 * 1024;
  static constexpr int STAGES_OFF = MT_HDR;
  static constexpr int TB = MT_BLOCKS * R * MC * 4;        // one fold buffer: [block][R][MC]
  static constexpr int TB_OFF = STAGES_OFF + NS * STAGE;
  static constexpr int BYTES = TB_OFF + 2 * TB;
  static constexpr int SMEM = BYTES + 1024;                // slack to align the base
  // the fold: each of the 32*TW fold threads owns FC columns of FRW rows
  static constexpr int FPT = R * MC / (32 * TW);           // (row, column) pairs per fold thread
  static constexpr int FC = FPT < MC ? FPT : MC;           // columns per fold thread
  static constexpr int FRW = FPT / FC;                     // rows per fold thread
  static constexpr int TPG = 32 * TW / (MC / FC);          // fold threads per column group
};

struct MtPlan {
  int tiles;     // row tiles x column chunks
  int CC;        // column chunks (of MC columns)
  int NSEG;      // segments per row (ceil(K / 512))
  const unsigned char* tabs;   // table records [CC][NSEG] in the workspace
};

// mbarriers in the header: stage full/empty, fold buffer full/empty
struct MtBars {
  uint64_t full[MT_NSMAX], empty[MT_NSMAX];
  uint64_t bfull[2], bempty[2];
};

// Untiled bulk copy global -> shared (16-byte aligned ends, a multiple of 16
// bytes), completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   sa(dst)),
               "l"(src), "r"(bytes), "r"(sa(bar))
               : "memory");
}

// The table of segment blockIdx.x for the column chunk blockIdx.y: the M = 1
// pipeline's scaled fp32 pairs of each column, side by side, and (fast mode)
// the block sums, in the record layout above.  Activations past M or K read
// as zero.  Exact form: step k of an item holds (code k of block 0, code k of
// block 1) * 2^-o(k); folded form: step 16*blk + CPW*p + j holds (code j of
// word 2p, of word 2p + 1) * 2^(FOLD_E - o(j)).  The block sums add the
// block's activations in the order of the dots (even and odd words serially,
// then together) and scale by 2^(b-1).
template <int BITS, bool FOLD, int MC, bool FUSED>
__global__ void __launch_bounds__(MT_TB_THREADS * MC)
    mt_table_kernel(const __half* x, const __half* r, const __half* gamma, float eps, __half* h_out, int M, int K,
                    int NSEG, unsigned char* tabs) {
  using RC = MtRec<MC>;
  constexpr int CPW = 32 / BITS, HALF = CPW / 2;
  __shared__ __align__(16) __half xs[2 * MC * 256];       // [half][m][256]
  __shared__ __align__(16) u64 rec[RC::TBLK / 8];
  extern __shared__ float nrm[];                           // fused: [MC][K/32] block sums, then [MC] inv
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // x (and r) come from the previous kernel, and it may still read the
  // workspace or h_out
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int s = blockIdx.x, m0 = blockIdx.y * MC, tt = threadIdx.x;
  for (int i = tt; i < RC::TBLK / 8; i += MT_TB_THREADS * MC) rec[i] = 0ull;
  if (FUSED) {
    // the residual add + RMSNorm of the fused definition, per column: warp
    // w takes column m0 + w, its lanes the block sums of squares of h =
    // fp16(x + r) (each serial over its 32 elements), lane 0 their serial
    // sum and inv = 1/sqrt(ss/K + eps) -- the same steps and order as the
    // M = 1 prologue, so the normalised activations are the same values
    const int NB = K / 32, w = tt >> 5, lane = tt & 31;
    float* bsum = nrm + w * NB;
    float* inv = nrm + MC * NB;
    if (m0 + w < M) {
      const __half* xc = x + (int64_t)(m0 + w) * K;
      const __half* rc = r + (int64_t)(m0 + w) * K;
      for (int b = lane; b < NB; b += 32) bsum[b] = block_sumsq(xc, rc, 32 * b, nullptr);
      __syncwarp();
      if (lane == 0) {
        float ss = 0.0f;
        for (int b = 0; b < NB; ++b) ss = __fadd_rn(ss, bsum[b]);
        inv[w] = rms_inv(ss, K, eps);
      }
    }
    __syncthreads();
  }
  for (int i = tt; i < MC * MT_KS / 8; i += MT_TB_THREADS * MC) {
    const int m = i / (MT_KS / 8), k = 8 * (i % (MT_KS / 8)), kk = s * MT_KS + k;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (m0 + m < M && kk < K) {
      const int64_t o = (int64_t)(m0 + m) * K + kk;
      if (FUSED) {
        // y = fp16((h * inv) * gamma), and h itself to h_out (this segment
        // of this chunk's columns)
        const uint4 xv = ldg16(reinterpret_cast<const uint4*>(x + o));
        const uint4 rv = ldg16(reinterpret_cast<const uint4*>(r + o));
        const uint4 gv = ldg16(reinterpret_cast<const uint4*>(gamma + kk));
        const float iv = nrm[MC * (K / 32) + m];
        uint16_t hh[8], yy[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const __half h = add_h(h_of(xv, e), h_of(rv, e));
          hh[e] = __half_as_ushort(h);
          yy[e] = __half_as_ushort(norm_h(h, iv, h_of(gv, e)));
        }
        memcpy(&v, yy, 16);
        if (h_out) {
          uint4 hv;
          memcpy(&hv, hh, 16);
          *reinterpret_cast<uint4*>(h_out + o) = hv;
        }
      } else {
        v = *reinterpret_cast<const uint4*>(x + o);
      }
    }
    *reinterpret_cast<uint4*>(xs + (k >> 8) * (MC * 256) + m * 256 + (k & 255)) = v;
  }
  __syncthreads();
  const int items = min(MT_ITEMS, (K - s * MT_KS) / 64);
  // 8 fp16 activations of column m from element k (a multiple of 8)
  auto chunk = [&](int m, int k, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(xs + (k >> 8) * (MC * 256) + m * 256 + (k & 255));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 h2 = u32_as_h2(w[e]);
      f[2 * e] = __low2float(h2);
      f[2 * e + 1] = __high2float(h2);
    }
  };
  // task (m, item, quarter): 8 steps of one item for one column, from two
  // 16-byte chunks of activations
  for (int task = tt; task < MC * items * 4; task += MT_TB_THREADS * MC) {
    const int m = task / (items * 4), iq = task % (items * 4), item = iq >> 2, q = iq & 3;
    const int hq = q & 1, blk = q >> 1;
    float A[8], Bv[8];
    if (!FOLD) {
      chunk(m, 64 * item + 8 * q, A);          // block 0, codes 8q ..
      chunk(m, 64 * item + 32 + 8 * q, Bv);    // block 1, codes 8q ..
    } else {
      const int a0 = 64 * item + 32 * blk + (BITS == 2 ? 8 : 16) * hq;
      chunk(m, a0, A);
      chunk(m, a0 + (BITS == 2 ? 16 : 8), Bv);
    }
    u64* dst = rec + (size_t)item * RC::TITEM + q * RC::OCT + m;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float v0, v1, sc;
      if (!FOLD) {
        sc = pow2f(-BITS * (((8 * q + i) % CPW) % HALF));
        v0 = A[i];
        v1 = Bv[i];
      } else {
        const int j = (8 * hq + i) % CPW;
        sc = pow2f(FOLD_E - BITS * (j % HALF));
        if (BITS == 8) {
          v0 = (i < 4) ? A[i] : Bv[i - 4];
          v1 = (i < 4) ? A[i + 4] : Bv[i];
        } else {
          v0 = A[i];
          v1 = Bv[i];
        }
      }
      dst[i * MC] = pk(__fmul_rn(v0, sc), __fmul_rn(v1, sc));
    }
  }
  if (FOLD) {
    float* ysum = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(rec) + RC::TAB);
    for (int task = tt; task < MC * 2 * items; task += MT_TB_THREADS * MC) {
      const int m = task / (2 * items), bl = task % (2 * items);
      float y[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float f[8];
        chunk(m, 32 * bl + 8 * c, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[8 * c + e] = f[e];
      }
      float S0 = 0.0f, S1 = 0.0f;
#pragma unroll
      for (int t16 = 0; t16 < 16; ++t16) {
        const int k0 = 2 * CPW * (t16 / CPW) + t16 % CPW;
        S0 = __fadd_rn(S0, y[k0]);
        S1 = __fadd_rn(S1, y[k0 + CPW]);
      }
      ysum[bl * MC + m] = __fmul_rn(__fadd_rn(S0, S1), (float)(1 << (BITS - 1)));
    }
  }
  __syncthreads();
  uint4* out = reinterpret_cast<uint4*>(tabs + ((size_t)blockIdx.y * NSEG + s) * RC::TBLK);
  for (int i = tt; i < RC::TBLK / 16; i += MT_TB_THREADS * MC) out[i] = reinterpret_cast<const uint4*>(rec)[i];
}

template <int BITS, bool FOLD, int U, int MC_>
__global__ void __launch_bounds__(MtLayout<BITS, U, MC_>::THREADS, 1)
    gemm_mt_kernel(GemvArgs a, MtPlan P, const __grid_constant__ CUtensorMap tm_codes,
                   const __grid_constant__ CUtensorMap tm_scales) {
  using L = MtLayout<BITS, U, MC_>;
  using RC = MtRec<MC_>;
  constexpr int R = L::R, MC = L::MC, CW = L::CW, UW = L::UW, NS = L::NS;
  constexpr int CPW = 32 / BITS, HALF = CPW / 2, WPB = 32 / CPW, NP = 16 / CPW;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  constexpr int CPI = BITS / 2;          // 16-byte chunks per item and row
  constexpr int IPB = 8 / CPI;           // items per 128-byte box
  static_assert((MC == 4 || MC == 8) && (L::FC == 8 || L::FC == 4 || L::FC == 2 || L::FC == 1) &&
                    R * MC == 32 * L::TW * L::FC * L::FRW && L::TPG * L::FRW == R,
                "tile shape");

  extern __shared__ unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((1024u - (sa(sm_raw) & 1023u)) & 1023u);
  MtBars* B = reinterpret_cast<MtBars*>(sm);
  volatile int* abort_f = reinterpret_cast<volatile int*>(sm + 512);
  int* err = &g_mt_error;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t perrow = a.perrow;

  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&B->full[s], 1);
      mbar_init(&B->empty[s], CW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B->bfull[b], CW);
      mbar_init(&B->bempty[b], L::TW);
    }
    *abort_f = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // the tables come from the table kernel, and the previous kernel may still
  // read y
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ------------------------------------------------------------ copies --
  if (warp == CW + L::TW) {
    if (lane == 0) {
      const uint32_t tx = (uint32_t)(L::NBOX * L::BOX + (perrow ? 0 : R * 32) + RC::TBLK);
      int g = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < P.tiles && !stop; t += gridDim.x) {
        const int r0 = (t / P.CC) * R, c = t % P.CC;
        const unsigned char* trec = P.tabs + (size_t)c * P.NSEG * RC::TBLK;
        for (int s = 0; s < P.NSEG; ++s, ++g) {
          const int slot = g % NS;
          if (g >= NS &&
              !mbar_wait_fast(&B->empty[slot], ((g / NS) - 1) & 1, abort_f, ERR_MT_TIMEOUT, err)) {
            stop = true;
            break;
          }
          if (*abort_f) {
            stop = true;
            break;
          }
          unsigned char* st = sm + L::STAGES_OFF + slot * L::STAGE;
          mbar_arrive_tx(&B->full[slot], tx);
#pragma unroll
          for (int b = 0; b < L::NBOX; ++b) tma_2d(st + b * L::BOX, &tm_codes, s * 8 * BITS + 16 * b, r0, &B->full[slot]);
          if (!perrow) tma_2d(st + L::SC_OFF, &tm_scales, s * 16, r0, &B->full[slot]);
          bulk_g2s(st + L::TBL_OFF, trec + (size_t)s * RC::TBLK, RC::TBLK, &B->full[slot]);
        }
      }
      // let every copy issued land before the CTA can exit
      for (int j = (g > NS ? g - NS : 0); j < g; ++j) mbar_drain(&B->full[j % NS], (j / NS) & 1, err);
    }
    return;
  }

  // --------------------------------------------------------- fold warps --
  if (warp >= CW) {
    // Thread tt owns FC columns of FRW rows of the tile (rows ri + TPG*k) and
    // adds each segment's block results in block order; after a tile's last
    // segment it stores the tile.
    constexpr int FC = L::FC, FRW = L::FRW, TPG = L::TPG;
    const int tt = tid - 32 * CW;   // 0 .. 32*L::TW - 1
    const int ri = tt % TPG, fc0 = (tt / TPG) * FC;
    float acc[FRW][FC];
#pragma unroll
    for (int k = 0; k < FRW; ++k)
#pragma unroll
      for (int c = 0; c < FC; ++c) acc[k][c] = 0.0f;
    int g = 0;
    for (int t = blockIdx.x; t < P.tiles; t += gridDim.x) {
      const int r0 = (t / P.CC) * R, m0 = (t % P.CC) * MC;
      for (int s = 0; s < P.NSEG; ++s, ++g) {
        const int bb = g & 1;
        const int items = min(MT_ITEMS, (a.K - s * MT_KS) / 64);
        if (!mbar_wait_fast(&B->bfull[bb], (g >> 1) & 1, abort_f, ERR_MT_TIMEOUT, err)) return;
#pragma unroll
        for (int k = 0; k < FRW; ++k) {
          const float* tb = reinterpret_cast<const float*>(sm + L::TB_OFF + bb * L::TB) + (ri + TPG * k) * MC + fc0;
#pragma unroll
          for (int bl = 0; bl < MT_BLOCKS; ++bl)
            if (bl < 2 * items) {
              if constexpr (FC == 8) {
                const float4 f = *reinterpret_cast<const float4*>(tb + bl * R * MC);
                const float4 f2 = *reinterpret_cast<const float4*>(tb + bl * R * MC + 4);
                acc[k][0] = __fadd_rn(acc[k][0], f.x);
                acc[k][1] = __fadd_rn(acc[k][1], f.y);
                acc[k][2] = __fadd_rn(acc[k][2], f.z);
                acc[k][3] = __fadd_rn(acc[k][3], f.w);
                acc[k][4] = __fadd_rn(acc[k][4], f2.x);
                acc[k][5] = __fadd_rn(acc[k][5], f2.y);
                acc[k][6] = __fadd_rn(acc[k][6], f2.z);
                acc[k][7] = __fadd_rn(acc[k][7], f2.w);
              } else if constexpr (FC == 4) {
                const float4 f = *reinterpret_cast<const float4*>(tb + bl * R * MC);
                acc[k][0] = __fadd_rn(acc[k][0], f.x);
                acc[k][1] = __fadd_rn(acc[k][1], f.y);
                acc[k][2] = __fadd_rn(acc[k][2], f.z);
                acc[k][3] = __fadd_rn(acc[k][3], f.w);
              } else if constexpr (FC == 2) {
                const float2 f = *reinterpret_cast<const float2*>(tb + bl * R * MC);
                acc[k][0] = __fadd_rn(acc[k][0], f.x);
                acc[k][1] = __fadd_rn(acc[k][1], f.y);
              } else {
                acc[k][0] = __fadd_rn(acc[k][0], tb[bl * R * MC]);
              }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B->bempty[bb]);
        if (s == P.NSEG - 1) {
#pragma unroll
          for (int k = 0; k < FRW; ++k) {
            const int64_t n = (int64_t)r0 + ri + TPG * k;
#pragma unroll
            for (int c = 0; c < FC; ++c) {
              const int col = m0 + fc0 + c;
              if (n < a.N && col < a.M) {
                float out = acc[k][c];
                if (perrow) out = __fadd_rn(0.0f, __fmul_rn(out, __half2float(a.scales[n])));
                const int64_t o = (int64_t)col * a.N + n;
                if (a.y_f16)
                  reinterpret_cast<__half*>(a.y)[o] = __float2half_rn(out);
                else
                  reinterpret_cast<float*>(a.y)[o] = out;
              }
              acc[k][c] = 0.0f;
            }
          }
        }
      }
    }
    return;
  }

  // ----------------------------------------------------- compute warps --
  bool ok = true;
  int g = 0;
  for (int t = blockIdx.x; t < P.tiles; t += gridDim.x) {
    for (int s = 0; s < P.NSEG; ++s, ++g) {
      const int slot = g % NS, b = g & 1;
      const int items = min(MT_ITEMS, (a.K - s * MT_KS) / 64);
      if (ok) ok = mbar_wait_fast(&B->full[slot], (g / NS) & 1, abort_f, ERR_MT_TIMEOUT, err);
      if (ok && g >= 2) ok = mbar_wait_fast(&B->bempty[b], ((g >> 1) - 1) & 1, abort_f, ERR_MT_TIMEOUT, err);

      // item `warp / CWI` of the segment for rows half `warp % CWI` of the
      // tile (lane: rows lane + 32 * (half * UW + u))
      const int item = warp / L::CWI, rh = (warp % L::CWI) * UW;
      if (ok && item < items) {
        const unsigned char* st = sm + L::STAGES_OFF + slot * L::STAGE;
        const u64* tabi = reinterpret_cast<const u64*>(st + L::TBL_OFF) + (size_t)item * RC::TITEM;
        const float* ysum = reinterpret_cast<const float*>(st + L::TBL_OFF + RC::TAB);
        float* tb = reinterpret_cast<float*>(sm + L::TB_OFF + b * L::TB);
        const unsigned char* cbox = st + (item / IPB) * L::BOX;
        const int ch0 = (item % IPB) * CPI;
        u64 wp[UW][BITS];   // the item's words as 64-bit pairs (2q, 2q + 1)
        uint32_t scw[UW];
#pragma unroll
        for (int u = 0; u < UW; ++u) {
          const int r = lane + 32 * (rh + u);
#pragma unroll
          for (int c = 0; c < CPI; ++c) {
            // 128-byte swizzle: chunk c of row r sits at chunk c ^ (r % 8)
            const ulonglong2 v =
                *reinterpret_cast<const ulonglong2*>(cbox + r * 128 + (((ch0 + c) ^ (lane & 7)) << 4));
            wp[u][2 * c] = v.x;
            wp[u][2 * c + 1] = v.y;
          }
          scw[u] = perrow ? 0u : *reinterpret_cast<const uint32_t*>(st + L::SC_OFF + r * 32 + item * 4);
        }
        if (FOLD) {
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            u64 acc2[UW][MC];
#pragma unroll
            for (int u = 0; u < UW; ++u)
#pragma unroll
              for (int mm = 0; mm < MC; ++mm) acc2[u][mm] = 0ull;
#pragma unroll
            for (int p = 0; p < NP; ++p) {
              u64 lo[UW], hi[UW];
#pragma unroll
              for (int u = 0; u < UW; ++u) {
                lo[u] = wp[u][blk * NP + p];
                hi[u] = lo[u] >> 16;
              }
#pragma unroll
              for (int j = 0; j < CPW; ++j) {
                const uint32_t m32 = MASK << (BITS * (j % HALF));
                const u64 mm64 = ((u64)m32 << 32) | m32;
                u64 v[UW];
#pragma unroll
                for (int u = 0; u < UW; ++u) v[u] = ((j < HALF) ? lo[u] : hi[u]) & mm64;
                const int tq = CPW * p + j;   // step 16*blk + tq
                const u64* yk = tabi + (2 * blk + (tq >> 3)) * RC::OCT + (tq & 7) * MC;
#pragma unroll
                for (int mm = 0; mm < MC; mm += 2) {
                  const ulonglong2 y2 = *reinterpret_cast<const ulonglong2*>(yk + mm);
#pragma unroll
                  for (int u = 0; u < UW; ++u) {
                    acc2[u][mm] = ffma2(y2.x, v[u], acc2[u][mm]);
                    acc2[u][mm + 1] = ffma2(y2.y, v[u], acc2[u][mm + 1]);
                  }
                }
              }
            }
            const int bl = 2 * item + blk;
            float bs[MC];
#pragma unroll
            for (int c4 = 0; c4 < MC; c4 += 4) {
              const float4 bS = *reinterpret_cast<const float4*>(ysum + bl * MC + c4);
              bs[c4] = bS.x;
              bs[c4 + 1] = bS.y;
              bs[c4 + 2] = bS.z;
              bs[c4 + 3] = bS.w;
            }
#pragma unroll
            for (int u = 0; u < UW; ++u) {
              const float sc = __half2float(__ushort_as_half((uint16_t)(blk ? (scw[u] >> 16) : (scw[u] & 0xFFFFu))));
              float o[MC];
#pragma unroll
              for (int mm = 0; mm < MC; ++mm) {
                float pe, po;
                upk(acc2[u][mm], pe, po);
                float pb = fold_block(__fadd_rn(pe, po), bs[mm]);
                if (!perrow) pb = __fmul_rn(pb, sc);
                o[mm] = pb;
              }
#pragma unroll
              for (int c4 = 0; c4 < MC; c4 += 4)
                *reinterpret_cast<float4*>(tb + (bl * R + lane + 32 * (rh + u)) * MC + c4) =
                    make_float4(o[c4], o[c4 + 1], o[c4 + 2], o[c4 + 3]);
            }
          }
        } else {
          uint32_t w[UW][2 * WPB];
#pragma unroll
          for (int u = 0; u < UW; ++u)
#pragma unroll
            for (int q = 0; q < BITS; ++q) {
              w[u][2 * q] = (uint32_t)wp[u][q];
              w[u][2 * q + 1] = (uint32_t)(wp[u][q] >> 32);
            }
          u64 acc2[UW][MC];
#pragma unroll
          for (int u = 0; u < UW; ++u)
#pragma unroll
            for (int mm = 0; mm < MC; ++mm) acc2[u][mm] = 0ull;
#pragma unroll
          for (int wi = 0; wi < WPB; ++wi) {
            uint32_t h0[UW], h1[UW];
#pragma unroll
            for (int u = 0; u < UW; ++u) {
              h0[u] = w[u][wi] >> 16;
              h1[u] = w[u][WPB + wi] >> 16;
            }
#pragma unroll
            for (int j = 0; j < CPW; ++j) {
              const int o = BITS * (j % HALF);
              const float offf = pow2f(23) + (float)(1 << (BITS - 1 + o));
              u64 v[UW];
#pragma unroll
              for (int u = 0; u < UW; ++u) {
                const uint32_t wa = (j < HALF) ? w[u][wi] : h0[u];
                const uint32_t wb = (j < HALF) ? w[u][WPB + wi] : h1[u];
                v[u] = decode2(wa, wb, MASK << o, pk(offf, offf));
              }
              const int tk = wi * CPW + j;   // step
              const u64* yk = tabi + (tk >> 3) * RC::OCT + (tk & 7) * MC;
#pragma unroll
              for (int mm = 0; mm < MC; mm += 2) {
                const ulonglong2 y2 = *reinterpret_cast<const ulonglong2*>(yk + mm);
#pragma unroll
                for (int u = 0; u < UW; ++u) {
                  acc2[u][mm] = ffma2(y2.x, v[u], acc2[u][mm]);
                  acc2[u][mm + 1] = ffma2(y2.y, v[u], acc2[u][mm + 1]);
                }
              }
            }
          }
#pragma unroll
          for (int u = 0; u < UW; ++u) {
            const float s_lo = __half2float(__ushort_as_half((uint16_t)(scw[u] & 0xFFFFu)));
            const float s_hi = __half2float(__ushort_as_half((uint16_t)(scw[u] >> 16)));
            const int r = lane + 32 * (rh + u);
            float o0[MC], o1[MC];
#pragma unroll
            for (int mm = 0; mm < MC; ++mm) {
              float p0, p1;
              upk(acc2[u][mm], p0, p1);
              o0[mm] = perrow ? p0 : __fmul_rn(p0, s_lo);
              o1[mm] = perrow ? p1 : __fmul_rn(p1, s_hi);
            }
#pragma unroll
            for (int c4 = 0; c4 < MC; c4 += 4) {
              *reinterpret_cast<float4*>(tb + ((2 * item) * R + r) * MC + c4) =
                  make_float4(o0[c4], o0[c4 + 1], o0[c4 + 2], o0[c4 + 3]);
              *reinterpret_cast<float4*>(tb + ((2 * item + 1) * R + r) * MC + c4) =
                  make_float4(o1[c4], o1[c4 + 1], o1[c4 + 2], o1[c4 + 3]);
            }
          }
        }
      }
      // the stage and this warp's share of the fold buffer are done
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&B->empty[slot]);
        mbar_arrive(&B->bfull[b]);
      }
    }
  }
}

}  // namespace

// ------------------------------------------------------------- launcher --

int read_mt_error(int clear, int* out) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_mt_error, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  if (clear && v) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_mt_error, &z, sizeof(int));
    if (e != cudaSuccess) return (int)e;
  }
  *out = v;
  return 0;
}

namespace {

// Launch on s, as a programmatic dependent of the previous kernel when PDL is
// on (every kernel here waits for its predecessor with griddepcontrol.wait).
template <typename... KArgs, typename... Args>
cudaError_t mt_launch(void (*kern)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t s,
                      Args... args) {
  if (pdl_enabled()) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
  }
  kern<<<grid, threads, smem, s>>>(args...);
  return cudaGetLastError();
}

size_t mt_table_bytes(int M, int K, int MC) {
  const size_t CC = (size_t)(M + MC - 1) / MC, NSEG = (size_t)(K + MT_KS - 1) / MT_KS;
  return CC * NSEG * (size_t)(MC == 8 ? MtRec<8>::TBLK : MtRec<4>::TBLK);
}

// The table kernel, then the tiles on its records (a.ws: the records).
template <int BITS, bool FOLD, int U, int MC>
int run_mt(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  using L = MtLayout<BITS, U, MC>;
  constexpr int R = L::R;
  auto kern = gemm_mt_kernel<BITS, FOLD, U, MC>;
  static thread_local KernCache cache;
  const DevInfo& d = dev_info();
  if ((size_t)L::SMEM > (size_t)d.max_smem_optin) return QMV_ERR_UNSUPPORTED;
  if (!a.ws || a.ws_bytes < mt_table_bytes(a.M, a.K, MC)) return QMV_ERR_WORKSPACE;
  int occ = 0;
  cudaError_t e = prep_kernel(kern, cache, L::THREADS, L::SMEM, &occ);
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  if (occ < 1) return QMV_ERR_UNSUPPORTED;
  // codes as UINT64 [N][row_bytes/8] (box 16 x R, 128-byte swizzle), scales
  // as UINT16 [N][K/32] (box 16 x R); rows past N are zero-filled
  const uint64_t row_bytes = (uint64_t)a.K * BITS / 8;
  CUtensorMap tmc, tms;
  if (!enc2d(&tmc, CU_TENSOR_MAP_DATA_TYPE_UINT64, a.codes, row_bytes / 8, (uint64_t)a.N, row_bytes, 16, R,
             CU_TENSOR_MAP_SWIZZLE_128B))
    return QMV_ERR_UNSUPPORTED;
  if (a.perrow)
    tms = tmc;   // unused
  else if (!enc2d(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.scales, (uint64_t)a.G, (uint64_t)a.N,
                  (uint64_t)a.G * 2, 16, R, CU_TENSOR_MAP_SWIZZLE_NONE))
    return QMV_ERR_UNSUPPORTED;
  MtPlan P;
  P.CC = (a.M + MC - 1) / MC;
  P.tiles = (int)(((int64_t)a.N + R - 1) / R) * P.CC;
  P.NSEG = (a.K + MT_KS - 1) / MT_KS;
  P.tabs = reinterpret_cast<const unsigned char*>(a.ws);
  if (a.fused) {
    // the fused residual add + RMSNorm runs in the table kernel
    const size_t nsm = ((size_t)MC * (a.K / 32) + MC) * sizeof(float);
    auto tk = mt_table_kernel<BITS, FOLD, MC, true>;
    if (nsm > 16 * 1024) e = cudaFuncSetAttribute(tk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)nsm);
    if (e == cudaSuccess)
      e = mt_launch(tk, dim3(P.NSEG, P.CC), MT_TB_THREADS * MC, nsm, s, a.x, a.r, a.gamma, a.eps, a.h_out, a.M, a.K,
                    P.NSEG, reinterpret_cast<unsigned char*>(a.ws));
  } else {
    e = mt_launch(mt_table_kernel<BITS, FOLD, MC, false>, dim3(P.NSEG, P.CC), MT_TB_THREADS * MC, 0, s, a.x,
                  (const __half*)nullptr, (const __half*)nullptr, 0.0f, (__half*)nullptr, a.M, a.K, P.NSEG,
                  reinterpret_cast<unsigned char*>(a.ws));
  }
  if (e == cudaSuccess) {
    const int grid = P.tiles < d.sms ? P.tiles : d.sms;
    e = mt_launch(kern, dim3(grid), L::THREADS, L::SMEM, s, a, P, tmc, tms);
  }
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  return QMV_OK;
}

// The tile shapes built: rows per lane U and columns MC.  8-column tiles
// share each code's mask between twice the paired FMAs; they fit shared
// memory with two ring stages, for int2 at U <= 4 and for int4 and int8 at
// U = 2.
struct MtChoice {
  int U, MC;
};
static bool mt_built(int bits, int U, int MC) {
  if (MC == 4) return U == 1 || U == 2 || (U == 4 && bits != 8);
  return U == 2 || (U == 4 && bits == 2);
}

// Estimated time of a tile shape, in SM cycles: whole rounds of tiles over
// the SMs, times the segments per tile, times the measured cost of one
// segment on GB300 (4 columns: about 4500 cycles for 128 rows, 2900 for 64,
// 32-row tiles priced on the same line; 8 columns: twice the paired FMAs at
// about 10 % better issue efficiency on the same fixed part).
static double mt_cost(int N, int M, int K, int U, int MC, int sms) {
  const int R = 32 * U;
  const int64_t tiles = (((int64_t)N + R - 1) / R) * ((M + MC - 1) / MC);
  const int64_t rounds = (tiles + sms - 1) / sms;
  const double seg = (MC == 4) ? 1300.0 + 25.0 * R : 1300.0 + 45.0 * R;
  return (double)rounds * ((K + MT_KS - 1) / MT_KS) * seg;
}

static MtChoice mt_choose(int N, int M, int K, int bits) {
  const int sms = dev_info().sms;
  MtChoice best{2, 4};
  double bc = mt_cost(N, M, K, 2, 4, sms);
  const MtChoice cand[] = {{4, 4}, {1, 4}, {2, 8}, {4, 8}};
  for (const MtChoice& c : cand) {
    if (!mt_built(bits, c.U, c.MC) || (c.MC == 8 && M < 5)) continue;
    const double t = mt_cost(N, M, K, c.U, c.MC, sms);
    if (t < bc) {
      bc = t;
      best = c;
    }
  }
  return best;
}

template <int BITS, bool FOLD>
int mt_bits(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  const MtChoice c = mt_choose(a.N, a.M, a.K, BITS);
  if (c.MC == 8) {
    if constexpr (BITS == 2)
      if (c.U == 4) return run_mt<BITS, FOLD, 4, 8>(a, s, err);
    return run_mt<BITS, FOLD, 2, 8>(a, s, err);
  }
  if (c.U == 1) return run_mt<BITS, FOLD, 1, 4>(a, s, err);
  if constexpr (BITS != 8)
    if (c.U == 4) return run_mt<BITS, FOLD, 4, 4>(a, s, err);
  return run_mt<BITS, FOLD, 2, 4>(a, s, err);
}

}  // namespace

static int launch_mtile_plain(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err);

size_t mt_workspace_bytes(int M, int N, int K, int bits, bool fused) {
  (void)fused;   // the fused residual add + RMSNorm needs no scratch of its own
  if (M < 2 || K % 256 != 0) return 0;
  const MtChoice c = mt_choose(N, M, K, bits);
  return mt_table_bytes(M, K, c.MC);
}

int launch_mtile(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err) {
  if (a.M < 2 || a.K % 256 != 0 || a.gather_rows || a.amax_ws) return QMV_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(a.x) & 15u) != 0) return QMV_ERR_UNSUPPORTED;
  if (!a.ws || a.ws_bytes < mt_workspace_bytes(a.M, a.N, a.K, bits, a.fused != 0)) return QMV_ERR_WORKSPACE;
  return launch_mtile_plain(a, bits, s, err);
}

static int launch_mtile_plain(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err) {
  if (a.folded) {
    switch (bits) {
      case 2: return mt_bits<2, true>(a, s, err);
      case 4: return mt_bits<4, true>(a, s, err);
      default: return mt_bits<8, true>(a, s, err);
    }
  }
  switch (bits) {
    case 2: return mt_bits<2, false>(a, s, err);
    case 4: return mt_bits<4, false>(a, s, err);
    default: return mt_bits<8, false>(a, s, err);
  }
}

}  // namespace qmv
