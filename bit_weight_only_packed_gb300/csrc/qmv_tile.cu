// qmv_tile.cu -- M-column tiles (2 <= M <= 32 token columns) on paired fp32
// arithmetic, for K a multiple of 64.
//
// What they compute ("raw-metal-loop-playbook", prefill-regimes table: keep
// each output scalar's K-dot in the single-token accumulation order and stage
// the weights across the M columns): every column of a tile is bit-identical
// to the M = 1 pipeline's result for that column, in both modes -- the exact
// form (the oracle's order) and the fast mode's folded-offset form (see
// qmv_decode.cuh), which the M = 1 pipeline also uses when K is a multiple of
// 256.
#include "qmv_prologue.cuh"

namespace qmv {

// ============================================ M-column tiles, paired fp32 ====
//
// The same computation as gemm_small_kernel for K a multiple of 64, on the
// arithmetic of the M = 1 pipeline: every 64-code item (two 32-code blocks)
// is decoded per position into the exact fp32 pair (v_k, v_{32+k}) * 2^o with
// two LOP3s and one paired subtract, and one fma.rn.f32x2 per column advances
// that column's two block chains, with the activations pre-scaled by 2^-o in
// shared memory ((y*2^-o)*(v*2^o) = y*v exactly, so each step is the oracle's
// rounded fp32 add).  With FOLD (fast mode) the masked fields are the
// operands, the activations are pre-scaled by 2^(FOLD_E - o) and each block
// is finished with its activation sum, as in the M = 1 pipeline.  Lanes are
// rows; warp w takes item w of each 512-code slab; a column's activation
// pairs are read as shared-memory broadcasts, two columns per 16-byte load;
// columns are processed 16 at a time.

constexpr int TL_WARPS = 8;
constexpr int TL_SLAB = TL_WARPS * 64;   // codes per slab
constexpr int TL_SB = TL_SLAB / 32;      // blocks per slab

template <int MT, int U> struct TileCfg {
  static constexpr int ROWS = 32 * U;                // rows per CTA (U per lane)
  static constexpr int PAIRS = ROWS * MT;
  static constexpr int PPT = (PAIRS + 255) / 256;
  static constexpr int MS = MT + 2;                  // padded column stride of the pair table
  static constexpr int YP = TL_WARPS * 32 * MS;      // activation pairs (u64) per slab
  static constexpr int TB = TL_SB * MT * ROWS;       // fold buffer floats
};

// Shared memory: activation pairs, fold buffer (also the fp16 staging of a
// slab), inv per column, the fused prologue's
// block sums of squares, and (FOLD) the slab's per-block activation sums.
template <int MT, int U>
__host__ __device__ inline size_t tile_smem_bytes(int NB, bool fused, bool fold) {
  using S = TileCfg<MT, U>;
  size_t b = (size_t)S::YP * 8 + (size_t)S::TB * 4 + (size_t)((MT + 3) & ~3) * 4;
  if (fused) b += (size_t)MT * NB * 4;
  if (fold) b += (size_t)MT * TL_SB * 4;
  return b;
}

template <int BITS, int MT, int U, bool FOLD>
__global__ void __launch_bounds__(256) gemm_tile_kernel(GemvArgs a) {
  using S = TileCfg<MT, U>;
  static_assert(MT % 2 == 0, "column chunks are whole pairs");
  constexpr int IW = 64 * BITS / 32;      // words per item
  constexpr int CPW = 32 / BITS, HALF = CPW / 2, WPB = 32 / CPW;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  constexpr int MTC = (MT < 16) ? MT : 16;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // blockIdx.y selects a chunk of MT token columns (column split when there
  // are few row tiles)
  const int mc0 = blockIdx.y * MT;
  a.x += (int64_t)mc0 * a.K;
  if (a.fused) {
    a.r += (int64_t)mc0 * a.K;
    if (a.h_out) a.h_out += (int64_t)mc0 * a.K;
  }
  a.y = a.y_f16 ? (void*)(reinterpret_cast<__half*>(a.y) + (int64_t)mc0 * a.N)
                : (void*)(reinterpret_cast<float*>(a.y) + (int64_t)mc0 * a.N);
  a.M = min(MT, a.M - mc0);
  const int K = a.K, NB = K / 32, M = a.M;
  const int64_t row0 = (int64_t)blockIdx.x * S::ROWS;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  u64* yp = reinterpret_cast<u64*>(smem_raw);                 // [item][k][m], stride MT+2
  float* tb = reinterpret_cast<float*>(yp + S::YP);           // [block][m][row]
  float* inv = tb + S::TB;
  float* bsum = inv + ((MT + 3) & ~3);
  float* ssl = bsum + (a.fused ? MT * NB : 0);   // FOLD: [m][TL_SB] 2^(b-1) * S

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

  for (int s0 = 0; s0 < K; s0 += TL_SLAB) {
    const int items = min(TL_WARPS, (K - s0) / 64);
    // stage the slab's activations: (1) coalesced 16-byte loads (the fused
    // path forms h and y here) into an fp16 buffer [m][512] that aliases the
    // fold buffer (free between the fold and the block sums); (2) re-layout
    // into fp32 pairs (y_k, y_{32+k}) * 2^-o(k), [item][k][m] with column
    // stride MT+2, threads walking k fastest (conflict-free reads and stores)
    __half* y16 = reinterpret_cast<__half*>(tb);
    for (int e = t; e < MT * items * 8; e += 256) {
      const int m = e / (items * 8), kk = 8 * (e % (items * 8));
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
      *reinterpret_cast<uint4*>(y16 + m * TL_SLAB + kk) = out;
    }
    __syncthreads();
    if (FOLD) {
      // block sums of the activations in the order of the dots (even and
      // odd words serially, then added), times 2^(b-1)
      for (int e = t; e < MT * 2 * items; e += 256) {
        const int m = e / (2 * items), bl = e % (2 * items);
        const __half* yb = y16 + m * TL_SLAB + 32 * bl;
        float S0 = 0.0f, S1 = 0.0f;
#pragma unroll
        for (int tt = 0; tt < 16; ++tt) {
          const int k0 = CPW * 2 * (tt / CPW) + tt % CPW;
          S0 = __fadd_rn(S0, __half2float(yb[k0]));
          S1 = __fadd_rn(S1, __half2float(yb[k0 + CPW]));
        }
        ssl[m * TL_SB + bl] = __fmul_rn(__fadd_rn(S0, S1), (float)(1 << (BITS - 1)));
      }
    }
    for (int e = t; e < items * 32 * MT; e += 256) {
      const int k = e & 31, m = (e >> 5) % MT, it = (e >> 5) / MT;
      const __half* yi = y16 + m * TL_SLAB + 64 * it;
      float v0, v1;
      if (!FOLD) {
        // step k: (code k of block 0, code k of block 1)
        const float sc = pow2f(-BITS * ((k % CPW) % HALF));
        v0 = __fmul_rn(__half2float(yi[k]), sc);
        v1 = __fmul_rn(__half2float(yi[32 + k]), sc);
      } else {
        // step k = 16*blk + CPW*p + j: (code j of word 2p, of word 2p + 1)
        const int blk = k >> 4, p = (k & 15) / CPW, j = (k & 15) % CPW;
        const float sc = pow2f(FOLD_E - BITS * (j % HALF));
        const int k0 = 32 * blk + CPW * 2 * p + j;
        v0 = __fmul_rn(__half2float(yi[k0]), sc);
        v1 = __fmul_rn(__half2float(yi[k0 + CPW]), sc);
      }
      yp[(it * 32 + k) * S::MS + m] = pk(v0, v1);
    }
    __syncthreads();

    if (FOLD && warp < items) {
      // folded form: item `warp` of this slab, one block at a time, for rows
      // lane + 32u of the tile; the words as 64-bit pairs (2q, 2q + 1)
      constexpr int NP = 16 / CPW;   // word pairs per block
      const int item = s0 / 64 + warp;
      u64 wp[U][IW / 2];
      uint32_t scw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t row = row0 + lane + 32 * u;
        scw[u] = 0u;
        if (row < a.N) {
          const ulonglong2* src =
              reinterpret_cast<const ulonglong2*>(a.codes + row * a.row_u4 + (int64_t)item * (IW / 4));
#pragma unroll
          for (int q = 0; q < IW / 4; ++q) {
            const ulonglong2 v = __ldg(src + q);
            wp[u][2 * q] = v.x;
            wp[u][2 * q + 1] = v.y;
          }
          if (!a.perrow) scw[u] = __ldg(reinterpret_cast<const unsigned int*>(a.scales + row * a.G + (int64_t)item * 2));
        } else {
#pragma unroll
          for (int q = 0; q < IW / 2; ++q) wp[u][q] = 0ull;
        }
      }
      const u64* yit = yp + (size_t)warp * 32 * S::MS;
#pragma unroll 1
      for (int c0 = 0; c0 < MT; c0 += MTC) {
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          u64 acc2[U][MTC];
#pragma unroll
          for (int u = 0; u < U; ++u)
#pragma unroll
            for (int mm = 0; mm < MTC; ++mm) acc2[u][mm] = 0ull;
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            u64 lo[U], hi[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              lo[u] = wp[u][blk * NP + p];
              hi[u] = lo[u] >> 16;
            }
#pragma unroll
            for (int j = 0; j < CPW; ++j) {
              const uint32_t m32 = MASK << (BITS * (j % HALF));
              const u64 mm64 = ((u64)m32 << 32) | m32;
              u64 v[U];
#pragma unroll
              for (int u = 0; u < U; ++u) v[u] = ((j < HALF) ? lo[u] : hi[u]) & mm64;
              const u64* yk = yit + (16 * blk + CPW * p + j) * S::MS + c0;
#pragma unroll
              for (int mm = 0; mm < MTC; mm += 2) {
                const ulonglong2 y2 = *reinterpret_cast<const ulonglong2*>(yk + mm);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                  acc2[u][mm] = ffma2(y2.x, v[u], acc2[u][mm]);
                  acc2[u][mm + 1] = ffma2(y2.y, v[u], acc2[u][mm + 1]);
                }
              }
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const float sc = __half2float(__ushort_as_half((uint16_t)(blk ? (scw[u] >> 16) : (scw[u] & 0xFFFFu))));
#pragma unroll
            for (int mm = 0; mm < MTC; ++mm) {
              float pe, po;
              upk(acc2[u][mm], pe, po);
              float pb = fold_block(__fadd_rn(pe, po), ssl[(c0 + mm) * TL_SB + 2 * warp + blk]);
              if (!a.perrow) pb = __fmul_rn(pb, sc);
              tb[((2 * warp + blk) * MT + c0 + mm) * S::ROWS + lane + 32 * u] = pb;
            }
          }
        }
      }
    } else if (!FOLD && warp < items) {
      // item `warp` of this slab for rows lane + 32u of the tile
      const int item = s0 / 64 + warp;
      uint32_t w[U][IW];
      float s_lo[U], s_hi[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t row = row0 + lane + 32 * u;
        uint32_t sc = 0u;
        if (row < a.N) {
          const uint4* src = a.codes + row * a.row_u4 + (int64_t)item * (IW / 4);
#pragma unroll
          for (int q = 0; q < IW / 4; ++q) {
            const uint4 v = ldg16(src + q);
            w[u][4 * q] = v.x; w[u][4 * q + 1] = v.y; w[u][4 * q + 2] = v.z; w[u][4 * q + 3] = v.w;
          }
          if (!a.perrow) sc = __ldg(reinterpret_cast<const unsigned int*>(a.scales + row * a.G + (int64_t)item * 2));
        } else {
#pragma unroll
          for (int q = 0; q < IW; ++q) w[u][q] = 0u;
        }
        s_lo[u] = __half2float(__ushort_as_half((uint16_t)(sc & 0xFFFFu)));
        s_hi[u] = __half2float(__ushort_as_half((uint16_t)(sc >> 16)));
      }
      const u64* yit = yp + (size_t)warp * 32 * S::MS;
#pragma unroll 1
      for (int c0 = 0; c0 < MT; c0 += MTC) {
        u64 acc2[U][MTC];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int mm = 0; mm < MTC; ++mm) acc2[u][mm] = 0ull;
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
            u64 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const uint32_t wa = (j < HALF) ? w[u][wi] : h0[u];
              const uint32_t wb = (j < HALF) ? w[u][WPB + wi] : h1[u];
              v[u] = decode2(wa, wb, MASK << o, pk(offf, offf));
            }
            const u64* yk = yit + (wi * CPW + j) * S::MS + c0;
#pragma unroll
            for (int mm = 0; mm < MTC; mm += 2) {
              const ulonglong2 y2 = *reinterpret_cast<const ulonglong2*>(yk + mm);
#pragma unroll
              for (int u = 0; u < U; ++u) {
                acc2[u][mm] = ffma2(y2.x, v[u], acc2[u][mm]);
                acc2[u][mm + 1] = ffma2(y2.y, v[u], acc2[u][mm + 1]);
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int mm = 0; mm < MTC; ++mm) {
            float p0, p1;
            upk(acc2[u][mm], p0, p1);
            const int r = lane + 32 * u;
            tb[((2 * warp) * MT + c0 + mm) * S::ROWS + r] = a.perrow ? p0 : __fmul_rn(p0, s_lo[u]);
            tb[((2 * warp + 1) * MT + c0 + mm) * S::ROWS + r] = a.perrow ? p1 : __fmul_rn(p1, s_hi[u]);
          }
      }
    }
    __syncthreads();

    // fold this slab's blocks, in order, into the (row, column) accumulators
    const int sbe = 2 * items;
#pragma unroll
    for (int i = 0; i < S::PPT; ++i) {
      const int pq = t + 256 * i;
      if (pq < S::PAIRS) {
        const int prow = pq % S::ROWS, pm = pq / S::ROWS;
        float v = acc[i];
        for (int b = 0; b < sbe; ++b) v = __fadd_rn(v, tb[(b * MT + pm) * S::ROWS + prow]);
        acc[i] = v;
      }
    }
    // the next slab's staging reuses the fold buffer
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < S::PPT; ++i) {
    const int pq = t + 256 * i;
    if (pq < S::PAIRS) {
      const int prow = pq % S::ROWS, pm = pq / S::ROWS;
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

// ============================================================ launcher ====

template <int BITS, int MT, int U>
static int run_tile(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  const int NB = a.K / 32;
  const bool fold = a.folded != 0;
  const size_t smem = tile_smem_bytes<MT, U>(NB, a.fused != 0, fold);
  const DevInfo& d = dev_info();
  if (smem > (size_t)d.max_smem_optin) return QMV_ERR_UNSUPPORTED;
  auto kern = fold ? gemm_tile_kernel<BITS, MT, U, true> : gemm_tile_kernel<BITS, MT, U, false>;
  static thread_local KernCache cache[2];
  cudaError_t e = prep_kernel(kern, cache[fold ? 1 : 0], 256, smem, nullptr);
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  const int64_t grid = ((int64_t)a.N + 32 * U - 1) / (32 * U);
  const int chunks = (a.M + MT - 1) / MT;
  kern<<<dim3((unsigned)grid, (unsigned)chunks), 256, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) { *err = e; return QMV_ERR_CUDA; }
  return QMV_OK;
}

// Two rows per lane (half the activation loads per FMA) where the registers
// and the fold buffer allow it; column chunk: the whole M, halved (down to 4)
// while there are fewer than 2 CTAs per SM of row tiles x chunks.
template <int BITS>
static int tile_bits(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  constexpr int U2 = (BITS == 8) ? 1 : 2;
  int mt = (a.M <= 4) ? 4 : (a.M <= 8) ? 8 : (a.M <= 16) ? 16 : 32;
  const int64_t sms2 = 2LL * dev_info().sms;
  while (mt > 4 && (((int64_t)a.N + 63) / 64) * ((a.M + mt - 1) / mt) < sms2) mt /= 2;
  if (mt == 4) return run_tile<BITS, 4, U2>(a, s, err);
  if (mt == 8) return run_tile<BITS, 8, U2>(a, s, err);
  if (mt == 16) return run_tile<BITS, 16, U2>(a, s, err);
  return run_tile<BITS, 32, 1>(a, s, err);
}

int launch_tile(const GemvArgs& a, int bits, cudaStream_t s, cudaError_t* err) {
  if (a.K % 64 != 0 || a.M < 1 || a.M > 32) return QMV_ERR_UNSUPPORTED;
  switch (bits) {
    case 2: return tile_bits<2>(a, s, err);
    case 4: return tile_bits<4>(a, s, err);
    default: return tile_bits<8>(a, s, err);
  }
}

}  // namespace qmv
