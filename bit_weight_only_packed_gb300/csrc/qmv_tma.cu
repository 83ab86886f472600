// qmv_tma.cu -- the M = 1 matvec as a warp-specialised pipeline (GB300).
//
// What it computes is exactly what the CUDA-core kernels compute (and the
// oracle): per output row, each 32-code block summed serially in k in fp32
// with exact products, scaled (group 32), and folded serially over blocks
// ("Gemma4 raw-Metal loop on A19", section "What moved the needle": int2 at
// 16 codes per word, exact products, fp32 in code order; the residual-add +
// RMSNorm fold into the matvec prologue).  Fast mode runs the folded-offset
// form of the same sums (qmv_decode.cuh).
//
// How (building blocks in qmv_pipe.cuh):
//   * Rows are processed in groups of R rows, each in NSEG segments of K.  A
//     producer warp moves each (group, segment) -- R rows of codes and their
//     group-32 scales -- into a ring of M1_NS shared-memory stages with two
//     2-D tensor copies completing on the stage's "full" mbarrier.  It runs
//     ahead of the math by up to M1_NS stages and starts before the prologue,
//     since weights do not depend on the activations.
//   * Compute warps: thread t owns one 64-code item (two 32-code blocks) of
//     RP rows in parallel, U rows after another, reading the item's
//     activations from a shared-memory table pre-scaled per bit offset.  Exact
//     form: a field becomes fp32 exactly by one LOP3 ((w & (mask << o)) |
//     0x4B000000 = 2^23 + u*2^o), one paired subtract gives v*2^o, and one
//     paired FMA advances both blocks' serial sums.  Folded form: one 64-bit
//     AND per field pair and one paired FMA.
//   * Block sums (scaled) go to a ring of M1_TB fold buffers; a dedicated
//     fold warp adds them serially per row (one lane per row) and writes y,
//     so the compute warps never wait at a CTA-wide barrier.
//   * Every mbarrier wait is bounded; on timeout the kernel records an error
//     code in the device error word, stops issuing, lets its own copies land
//     and returns.
#include "qmv_pipe.cuh"

namespace qmv {

__device__ int g_qmv_error = 0;

using namespace pipe;

// Copy-ring stages and fold buffers of this kernel: three of each (against
// four stages and two fold buffers: the decode layer 923.6 -> 934.8 GB/s and
// the int4 262144 x 5376 lm_head 4.82 -> 4.94 TB/s) -- a third fold buffer
// lets the compute warps run two stages ahead of the fold warp, and the
// smaller ring pays for it in shared memory.
constexpr int M1_NS = 3, M1_TB = 3;
static_assert(8 * (2 * M1_NS + 2 * M1_TB) <= 96, "the kernel's mbarriers end below its flags at byte 96");

template <int BITS, bool PERROW, bool FUSED, bool EXACT, int U, int MAXT>
__global__ void __launch_bounds__(MAXT, (MAXT <= 320) ? 2 : 1)
    gemv_tma_kernel(GemvArgs a, TmaPlan P, const __grid_constant__ CUtensorMap tm_codes,
                    const __grid_constant__ CUtensorMap tm_scales) {
  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);
  uint64_t* empty = full + M1_NS;
  uint64_t* tfull = empty + M1_NS;
  uint64_t* tempty = tfull + M1_TB;
  volatile int* abort_f = reinterpret_cast<volatile int*>(sm + 96);
  float* inv_sh = reinterpret_cast<float*>(sm + 100);
  float* y2f = reinterpret_cast<float*>(sm + P.y_off);     // activation table
  float* ysum = reinterpret_cast<float*>(sm + P.ysum_off); // folded form: 2^(b-1) * S per block
  unsigned char* stages = sm + P.stage_off;
  float* tbuf = reinterpret_cast<float*>(sm + P.tbuf_off);
  int* ids_sh = reinterpret_cast<int*>(sm + P.ids_off);   // expert gather: selected ids
  int* err = &g_qmv_error;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = P.R;
  const int GS = P.KS / 32 + 4;          // fold-buffer row stride (16-byte aligned rows)
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
    if (threadIdx.x == 0) atomicCAS(err, 0, ERR_SMEM_ALIGN);
    return;
  }
  if (threadIdx.x == 0) {
    // consumers arrive once per warp (lane 0, after __syncwarp orders the
    // lanes' shared-memory accesses before its release)
    for (int s = 0; s < M1_NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], P.Tc / 32);
    }
    for (int b = 0; b < M1_TB; ++b) {
      mbar_init(&tfull[b], P.Tc / 32);
      mbar_init(&tempty[b], 1);
    }
    *abort_f = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ------------------------------------------------------------ producer --
  if (warp == 0) {
    if (a.gather_rows) {
      // the expert ids may come from the previous kernel: wait for it, then
      // keep them in shared memory (the fold warp reads them there, after
      // the stage barriers that follow these stores)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int t = lane; t < a.gather_n; t += 32) ids_sh[t] = a.gather_ids[t];
      __syncwarp();
    }
    int issued = 0;
    int seg = 0;
    int64_t g = blockIdx.x;
    for (int i = 0; i < my_stages; ++i) {
      const int s = i % M1_NS;
      if (i >= M1_NS && !mbar_wait_fast(&empty[s], ((i / M1_NS) - 1) & 1, abort_f, ERR_TIMEOUT_EMPTY, err)) break;
      if (*abort_f) break;
      const int64_t r0 = group_rows(a, R, g, ids_sh).phys0;
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
      for (int j = (issued > M1_NS ? issued - M1_NS : 0); j < issued; ++j)
        mbar_drain(&full[j % M1_NS], (j / M1_NS) & 1, err);
    return;
  }

  // ------------------------------------------- prologue (warps 1 .. end) --
  // Activations, residual and gamma may come from the previous kernel, and
  // the outputs may still be read by it: wait for it to complete (no-op
  // without a programmatic launch).  The producer above never waits: packed
  // weights are not written by the kernels a matvec overlaps.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the fold buffer is free until the main loop: it holds the block sums
  build_table<BITS, FUSED, EXACT>(a, y2f, ysum, tbuf, inv_sh, (blockIdx.x == 0) ? a.h_out : nullptr,
                                  threadIdx.x - 32, 32 + P.Tc, 1);
  named_bar(1, 32 + P.Tc);

  // ---------------------------------------------------------- fold warp --
  if (warp == 1) {
    float acc = 0.0f;   // this lane's row: group-32 accumulator, or the per-row block sum
    unsigned long long best = 0ull;   // argmax epilogue: this lane's best key
    int seg = 0;
    int64_t g = blockIdx.x;
    for (int i = 0; i < my_stages; ++i) {
      const int tb = i % M1_TB;
      if (!mbar_wait_fast(&tfull[tb], (i / M1_TB) & 1, abort_f, ERR_TIMEOUT_TFULL, err)) break;
      const GroupRows gr = group_rows(a, R, g, ids_sh);
      if (!gr.ok && lane == 0 && seg == 0) atomicCAS(err, 0, ERR_BAD_EXPERT);
      fold_stage(a, P, tbuf + (size_t)tb * R * GS, GS, lane, gr, seg, acc, a.amax_ws ? &best : nullptr);
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[tb]);
      if (++seg == P.NSEG) {
        seg = 0;
        g += gridDim.x;
      }
    }
    if (a.amax_ws) amax_finish(a, best, lane);
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
    const int s = i % M1_NS;
    const int tb = i % M1_TB;
    if (!mbar_wait_fast(&full[s], (i / M1_NS) & 1, abort_f, ERR_TIMEOUT_FULL, err)) break;
    if (i >= M1_TB && !mbar_wait_fast(&tempty[tb], ((i / M1_TB) - 1) & 1, abort_f, ERR_TIMEOUT_TEMPTY, err)) break;
    const int rows = a.gather_rows ? group_rows(a, R, g, ids_sh).rows
                                   : (int)min((int64_t)R, (int64_t)a.N - g * R);
    if (active)
      compute_stage<BITS, PERROW, EXACT, U>(stages + (size_t)s * P.stage_bytes, P, c, rp, seg, rows, y2s,
                                            ysum, tbuf + (size_t)tb * R * GS, GS);
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

// Plan for about `tc_target` compute threads and U rows per thread
// (RP*U <= 32 rows per group: one fold lane per row), in segments of at most
// ks_max codes.
static bool tma_plan(int N, int K, int bits, bool perrow, int tc_target, int U, TmaPlan* P,
                     int ks_max = 2048) {
  if (K % 256 != 0) return false;
  const int KS = tma_segment(K, ks_max);
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
  P->tbuf_off = tma_round16(P->stage_off + M1_NS * P->stage_bytes);
  {
    const int fold = M1_TB * P->R * (P->KS / 32 + 4) * 4;
    const int bsum = (K / 32) * 4;
    P->ids_off = P->tbuf_off + tma_round16(fold > bsum ? fold : bsum);
  }
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
// (K_seg / 32) x R.  tensor_maps caches them per thread (a few entries).
bool encode_pack_maps(const GemvArgs& a, const TmaPlan& P, CUtensorMap* tc, CUtensorMap* ts) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)(P.row_bytes / 8), (cuuint64_t)a.N};
    const cuuint64_t strides[1] = {(cuuint64_t)P.row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(P.seg_bytes / 8), (cuuint32_t)P.R};
    const cuuint32_t es[2] = {1, 1};
    if (enc(tc, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, (void*)a.codes, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  if (a.perrow) {
    *ts = *tc;   // unused
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 32), (cuuint64_t)a.N};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 32) * 2};
    const cuuint32_t box[2] = {(cuuint32_t)(P.KS / 32), (cuuint32_t)P.R};
    const cuuint32_t es[2] = {1, 1};
    if (enc(ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (void*)a.scales, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

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
  Entry e;
  e.codes = a.codes;
  e.scales = a.scales;
  e.N = a.N;
  e.K = a.K;
  e.bits = bits;
  e.R = P.R;
  e.KS = P.KS;
  if (!encode_pack_maps(a, P, &e.c, &e.s)) return false;
  cache[next] = e;
  next = (next + 1) % 8;
  if (valid < 8) ++valid;
  *tc = e.c;
  *ts = e.s;
  return true;
}

// Shared memory of a plan: up to the fold buffer (2 x R rows x (KS/32 + 1)
// floats, which also holds the fused prologue's K/32 block sums before the
// main loop), then room for GATHER_MAX expert ids.
static size_t tma_smem(const TmaPlan& P, int /*K*/) {
  return (size_t)P.ids_off + (size_t)GATHER_MAX * 4;
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
    if (U == 2) return run_tma<BITS, PERROW, FUSED, EXACT, 2, 576>(a, P, s, err, occ_only);
    if (U == 1) return run_tma<BITS, PERROW, FUSED, EXACT, 1, 576>(a, P, s, err, occ_only);
    return QMV_ERR_UNSUPPORTED;
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
// least 3 row groups per CTA slot when N allows it (load balance).  A small
// matrix (fewer than two such groups per CTA slot) may instead take the
// ~512-thread plan with one row per thread, when that shortens the busiest
// slot (ceil(groups / slots) stages, each a fixed part plus R rows).  The
// choice is cached per shape.
template <int BITS>
static int tma_bits(const GemvArgs& a, cudaStream_t s, cudaError_t* err) {
  struct Key { int N, K, perrow, fused, folded, gather, dev; };
  struct Entry { Key k; TmaPlan p; bool ok; };
  static thread_local Entry cache[16];
  static thread_local int next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  // rows the launch covers: the pack's, or the selected experts' (gather)
  const int Nl = a.gather_rows ? a.gather_n * a.gather_rows : a.N;
  auto gather_groups = [&](TmaPlan P) {
    if (a.gather_rows) P.ngroups = a.gather_n * ((a.gather_rows + P.R - 1) / P.R);
    return P;
  };
  const Key key{Nl, a.K, a.perrow, a.fused, a.folded, a.gather_rows, dev};
  for (int i = 0; i < 16; ++i) {
    const Key& k = cache[i].k;
    if (cache[i].ok && k.N == key.N && k.K == key.K && k.perrow == key.perrow &&
        k.fused == key.fused && k.folded == key.folded && k.gather == key.gather && k.dev == key.dev)
      return tma_dispatch<BITS>(a, gather_groups(cache[i].p), s, err, nullptr);
  }
  const int sms = dev_info().sms;
  TmaPlan best{};
  int best_score = -1;
  // small matrices (fewer than two full groups per CTA slot): a plan with
  // half-size groups (16 rows) -- one row per thread on 512 compute threads,
  // or, when K spans six or more segments, two rows per thread on 256 --
  // spreads the rows over more CTAs; it is taken when its busiest slot has
  // less to do.  Measured under graphs with programmatic dependent launch:
  // two rows per thread amortise each of many stages better (down
  // 2048x16384 int2 in a 30-layer token: 977 against 928 tok/s for the
  // token), while with up to four segments the 512-thread CTA is faster
  // (down 2048x8192 int2 in the decode layer: 22.75 against 23.65 us)
  TmaPlan small{};
  int64_t small_cost = -1, best_slots = 1;
  for (int tc : {256, 512}) {
    for (int U : {4, 2, 1}) {
      if (BITS == 8 && U > 2) continue;
      if (tc > 256 && U > 2) continue;
      if (tc <= 256 && U < 2) continue;
      TmaPlan P;
      if (!tma_plan(Nl, a.K, BITS, a.perrow != 0, tc, U, &P)) continue;
      if (tma_smem(P, a.K) > (size_t)dev_info().max_smem_optin) continue;
      int occ = 0;
      if (tma_dispatch<BITS>(a, gather_groups(P), s, err, &occ) != QMV_OK || occ < 1) continue;
      const TmaPlan Pg = gather_groups(P);
      const int64_t slots = (int64_t)occ * sms;
      const int64_t cost = ((Pg.ngroups + slots - 1) / slots) * (16 + P.R);
      if (U == 1 || (U == 2 && tc == 256 && P.R <= 16 && P.NSEG >= 6)) {
        if (small_cost < 0 || cost < small_cost || (cost == small_cost && U == 2)) {
          small_cost = cost;
          small = P;
        }
        if (U == 1) continue;
      }
      int score = occ * (P.Tc / 32) * 64 + P.R;
      // int4 is bound by the activation-table loads, which four rows per lane
      // halve: on large int4 matrices that beats a second CTA per SM (one
      // CTA of 224 compute threads at U = 4 against two of 256 at U = 2 on
      // the 262144 x 5376 lm_head: 4.82 against 4.24 TB/s)
      if (BITS == 4 && U == 4) score += 16 * 64;
      if ((int64_t)Pg.ngroups < 3LL * occ * sms && U > 2) score -= 64 * 64;   // balance
      if (score > best_score) {
        best_score = score;
        best = P;
        best_slots = slots;
      }
    }
  }
  if (best_score < 0) return QMV_ERR_UNSUPPORTED;
  if (small_cost >= 0) {
    const TmaPlan Bg = gather_groups(best);
    const int64_t best_cost = ((Bg.ngroups + best_slots - 1) / best_slots) * (16 + best.R);
    if ((int64_t)Bg.ngroups < 2 * best_slots && small_cost < best_cost) best = small;
  }
  // few rows over a long K (at most one 16-row group per SM): segments of
  // 4096 codes and four rows per thread on 256 compute threads, which halves
  // the activation-table reads per code against two rows per thread.
  // Measured on the int2 down projection 2048 x 16384 of a 30-layer decode
  // token (graphs with programmatic dependent launch): 877.5 -> 858.9 us a
  // token; 16 compute warps at two rows per thread gain nothing.
  if (BITS != 8 && a.K >= 16384 && a.K % 4096 == 0) {
    TmaPlan P;
    int occ = 0;
    if (tma_plan(Nl, a.K, BITS, a.perrow != 0, 256, 4, &P, 4096) && P.R == 16 &&
        tma_smem(P, a.K) <= (size_t)dev_info().max_smem_optin &&
        tma_dispatch<BITS>(a, gather_groups(P), s, err, &occ) == QMV_OK && occ >= 1 &&
        (int64_t)gather_groups(P).ngroups <= (int64_t)sms)
      best = P;
  }
  cache[next] = Entry{key, best, true};
  next = (next + 1) % 16;
  return tma_dispatch<BITS>(a, gather_groups(best), s, err, nullptr);
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
int read_chain_error(int clear, int* out);
int read_mt_error(int clear, int* out);

int read_device_error(int clear, int* out) {
  int t = 0, ch = 0, mt = 0;
  const int et = read_tc_error(clear, &t);
  if (et != 0) return et;
  const int ec = read_chain_error(clear, &ch);
  if (ec != 0) return ec;
  const int em = read_mt_error(clear, &mt);
  if (em != 0) return em;
  if (mt) t = mt;
  if (ch) t = ch;
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
